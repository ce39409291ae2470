"""GPU test of tq_attn_decode_noalloc, the decode entry point for callers that cannot
allocate device memory at decode time (frozen memory pools, plugins whose host framework
forbids cudaMalloc during a request): it must give the same outputs as tq_attn_decode with
a caller-provided workspace, on two calls in a row (the static scratch keeps the previous
call's contents), and reject requests larger than its 4 MiB scratch.

The file name makes pytest collect it last."""
import ctypes

import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import binding

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("d,b,G", [(128, 3, 4), (128, 3, 16), (64, 2, 2)])
def test_noalloc_matches_workspace_decode(d, b, G):
    B, H, T = 2, 2, 700
    ctx = tq.Context(d, b, seed=3)
    cache = ctx.alloc_cache(B, H, T)
    gen = torch.Generator().manual_seed(11)
    k = torch.randn(B, H, T, d, generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, T, d, generator=gen).to(torch.bfloat16).cuda()
    ctx.quantize_kv(k, v, torch.zeros(B, dtype=torch.int32, device="cuda"), cache, T)
    lens = torch.tensor([T, 301], dtype=torch.int32, device="cuda")
    ws = ctx.alloc_workspace(B, G * H, H, T)
    for call in range(2):
        q = torch.randn(B, G * H, d, generator=gen).cuda()
        ref = torch.empty_like(q)
        ctx.attn_decode(q, cache, lens, H, T, ref, ws)
        got = torch.full_like(q, float("nan"))
        rc = binding.tq_attn_decode_noalloc(ctx.handle, _ptr(q), B, G * H, H, _ptr(cache), _ptr(lens), T, _ptr(got),
                                            None, _stream())
        assert rc == tq.TQ_OK, tq.tq_status_string(rc)
        assert ctx.device_status() == tq.TQ_OK
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.isfinite(g)), call
        # the same kernels on the same inputs: identical up to the parity bar of the suite
        assert np.linalg.norm(g - r) <= 1e-6 * np.linalg.norm(r), call
    ctx.close()


def test_noalloc_rejects_requests_beyond_its_scratch():
    ctx = tq.Context(128, 3, seed=0)
    need = ctx.workspace_bytes(64, 1024, 64, 1 << 20)
    assert need > (4 << 20)
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    lens = torch.zeros(64, dtype=torch.int32, device="cuda")
    rc = binding.tq_attn_decode_noalloc(ctx.handle, _ptr(dummy), 64, 1024, 64, _ptr(dummy), _ptr(lens), 1 << 20,
                                        _ptr(dummy), None, _stream())
    assert rc == tq.TQ_ESCRATCH
    ctx.close()


def test_noalloc_returns_the_same_errors_as_decode():
    """A call the forced kernel cannot serve (the e2m1 tcgen05 kernel takes at most 8 query
    heads per KV head; here 12) and a group size that does not divide give tq_attn_decode's own
    error codes, not a generic one."""
    B, H, T, d = 1, 2, 256, 128
    ctx = tq.Context(d, 3, seed=0)
    ctx.set_decode_path("tc4")
    cache = ctx.alloc_cache(B, H, T)
    q = torch.zeros(B, 24, d, device="cuda")
    out = torch.empty_like(q)
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    rc_ref = binding.tq_attn_decode(ctx.handle, _ptr(q), B, 24, H, _ptr(cache), _ptr(lens), T, _ptr(out), None,
                                    _ptr(ws), ws.numel(), _stream())
    rc = binding.tq_attn_decode_noalloc(ctx.handle, _ptr(q), B, 24, H, _ptr(cache), _ptr(lens), T, _ptr(out), None,
                                        _stream())
    assert rc == rc_ref == tq.TQ_EUNSUPPORTED
    q3 = torch.zeros(B, 6, d, device="cuda")          # 6 query heads over 4 KV heads
    rc = binding.tq_attn_decode_noalloc(ctx.handle, _ptr(q3), B, 6, 4, _ptr(cache), _ptr(lens), T, _ptr(q3), None,
                                        _stream())
    assert rc == tq.TQ_EINVAL
    ctx.close()
