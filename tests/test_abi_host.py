"""CPU checks of the C-ABI library: it loads, exports every declared entry point, its host
argument checks reject bad input without touching a GPU, and its host-side set-up (seeded
Pi and S, Lloyd-Max codebooks) matches the oracle's independent implementation."""
import ctypes

import numpy as np
import pytest

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import binding
from oracle import codebook as ocb
from oracle import rotation as orot


def test_library_exports_every_declared_function():
    names = binding.header_functions()
    assert len(names) >= 13
    L = tq.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert missing == []
    assert set(binding._SIGS) == set(names)


def test_status_strings():
    assert tq.tq_status_string(0) == "ok"
    for code in range(-8, 0):
        assert tq.tq_status_string(code) != "unknown status"


@pytest.mark.parametrize("d", [8, 64, 128, 256])
def test_rotation_matches_oracle(d):
    pi = np.array(tq.tq_make_rotation(d, 0)).reshape(d, d)
    ref = orot.haar_rotation(d, 0)
    assert np.max(np.abs(pi - ref)) <= 1e-12
    assert np.max(np.abs(pi.T @ pi - np.eye(d))) <= 1e-12


@pytest.mark.parametrize("seed", [0, 1, 12345])
def test_projection_matches_oracle(seed):
    s = np.array(tq.tq_make_projection(128, 128, seed)).reshape(128, 128)
    ref = orot.qjl_matrix(128, 128, seed)
    assert np.max(np.abs(s - ref)) <= 1e-12


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("levels", [2, 4, 8, 16, 32])
def test_codebook_matches_oracle(d, levels):
    c, t = tq.tq_make_codebook(d, levels)
    rc, rt = ocb.codebook(d, levels)
    assert np.max(np.abs(np.array(c) - rc)) <= 1e-12
    assert np.max(np.abs(np.array(t) - rt)) <= 1e-12
    assert t[levels // 2 - 1] == 0.0


def test_host_argument_checks_need_no_gpu():
    L = tq.lib()
    out = ctypes.c_void_p()
    assert L.tq_ctx_create(100, 3, 100, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_create(128, 6, 128, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_create(128, 3, 64, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_create(128, 3, 128, 0, 0, None) == tq.TQ_EINVAL
    assert L.tq_quantize_kv(None, None, None, 1, 1, 1, None, None, 1, None) == tq.TQ_EINVAL
    assert L.tq_attn_decode(None, None, 1, 1, 1, None, None, 1, None, None, None, 0, None) == tq.TQ_EINVAL
    assert L.tq_cache_bytes(None, 1, 1, 1) == 0
    assert L.tq_decode_workspace_bytes(None, 1, 1, 1, 1) == 0
    assert L.tq_get_device_status(None, None) == tq.TQ_EINVAL
    assert L.tq_ctx_set_decode_path(None, tq.TQ_DECODE_TC) == tq.TQ_EINVAL
    c = (ctypes.c_double * 4)()
    assert L.tq_make_codebook(2, 4, c, c) == tq.TQ_EINVAL
    assert L.tq_make_codebook(128, 65, c, c) == tq.TQ_EINVAL


def test_host_argument_checks_of_the_extension_calls():
    """Format version 2, Sparse V, strided input, the paged pool and the scan reject bad
    arguments on the host (no GPU needed)."""
    L = tq.lib()
    out = ctypes.c_void_p()
    # format version 2: widths 1..5, d in {64, 128, 256}
    assert L.tq_ctx_create_kv(128, 7, 3, 1, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_create_kv(128, 3, 0, 0, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_create_kv(96, 3, 3, 1, 0, 0, ctypes.byref(out)) == tq.TQ_EUNSUPPORTED
    assert L.tq_ctx_set_sparse_v(None, 0.1) == tq.TQ_EINVAL
    st = (ctypes.c_int64 * 6)(0, 0, 128, 0, 0, 128)
    assert L.tq_quantize_kv_strided(None, None, None, st, 1, 1, 1, None, None, 1, None) == tq.TQ_EINVAL
    assert L.tq_quantize_kv_strided(None, None, None, None, 1, 1, 1, None, None, 1, None) == tq.TQ_EINVAL
    # paged pool: a missing pool or table, no blocks or no table columns
    assert L.tq_paged_pool_bytes(None, 1, 1) == 0
    assert L.tq_quantize_kv_paged(None, None, None, 1, 1, 1, None, None, 1, None, 1, None) == tq.TQ_EINVAL
    assert L.tq_quantize_kv_paged_strided(None, None, None, st, 1, 1, 1, None, None, 1, None, 1, None) == tq.TQ_EINVAL
    assert L.tq_attn_decode_paged(None, None, 1, 1, 1, None, 1, None, 1, None, None, None, None, 0,
                                  None) == tq.TQ_EINVAL
    assert L.tq_dequantize_kv_paged(None, None, 1, None, 1, 1, 1, None, 1, None, None, None) == tq.TQ_EINVAL
    # scan
    assert L.tq_ip_topk_workspace_bytes(None, 1, 1, 1, 1) == 0
    assert L.tq_ip_topk(None, None, 1, 1, 1, None, None, 1, 10, None, None, None, 0, None) == tq.TQ_EINVAL
    assert L.tq_ip_topk_paged(None, None, 1, 1, 1, None, 1, None, 1, None, 10, None, None, None, 0,
                              None) == tq.TQ_EINVAL


def test_binding_reads_strides_of_a_token_major_view():
    import torch
    B, T, H, d = 2, 5, 3, 128
    k = torch.zeros(B, T, H, d, dtype=torch.bfloat16)
    view = k.permute(0, 2, 1, 3)   # the quantizer's [B, H, T, d] view of a projection output
    st = tq.Context._kv_strides(view, view)
    assert list(st) == [T * H * d, d, H * d] * 2
    with pytest.raises(tq.TQError):
        tq.Context._kv_strides(view.transpose(2, 3), view.transpose(2, 3))   # d not contiguous
