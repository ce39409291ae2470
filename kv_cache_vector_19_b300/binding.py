"""ctypes binding of ``libtq.so``: the same entry points as ``include/tq.h``.

Argument marshalling only.  Every step of the quantize / decode path runs in the library's
CUDA kernels; PyTorch is used here for nothing but device memory and the current stream.
If the shared library cannot be built or loaded, every call raises: there is no fallback.
"""
import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "tq.h")
LIB_PATH = os.path.join(PKG, "libtq.so")

TQ_OK = 0
TQ_EINVAL = -1
TQ_EUNSUPPORTED = -2
TQ_ECUDA = -3
TQ_ETIMEOUT = -4
TQ_EBOUNDS = -5
TQ_ENOMEM = -6
TQ_ENOTCONV = -7
TQ_ESCRATCH = -8
TQ_TOPK_MAX = 1024
TQ_DECODE_AUTO, TQ_DECODE_SIMT, TQ_DECODE_MMA, TQ_DECODE_TC, TQ_DECODE_TC4 = 0, 1, 2, 3, 4
DECODE_PATHS = {"auto": TQ_DECODE_AUTO, "simt": TQ_DECODE_SIMT, "mma": TQ_DECODE_MMA, "tc": TQ_DECODE_TC,
                "tc4": TQ_DECODE_TC4}
PAGE_TOKENS = 128
# kernels one call launches (the benchmark reports launch counts from these)
QUANTIZE_LAUNCHES = 1
DECODE_LAUNCHES = 3

_lock = threading.Lock()
_lib = None

_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_dp = ctypes.POINTER(ctypes.c_double)

# name -> (restype, argtypes)
_SIGS = {
    "tq_make_codebook": (_c_int, [_c_int, _c_int, _dp, _dp]),
    "tq_make_rotation": (_c_int, [_c_int, ctypes.c_uint64, _dp]),
    "tq_make_projection": (_c_int, [_c_int, _c_int, ctypes.c_uint64, _dp]),
    "tq_ctx_create": (_c_int, [_c_int, _c_int, _c_int, ctypes.c_uint64, _c_int, ctypes.POINTER(_vp)]),
    "tq_ctx_create_kv": (_c_int, [_c_int, _c_int, _c_int, _c_int, ctypes.c_uint64, _c_int, ctypes.POINTER(_vp)]),
    "tq_ctx_destroy": (None, [_vp]),
    "tq_page_bytes": (_c_size, [_vp]),
    "tq_cache_bytes": (_c_size, [_vp, _c_int, _c_int, _c_int]),
    "tq_ctx_get_constants": (_c_int, [_vp, _dp, _dp, _dp, _dp, _dp, _dp]),
    "tq_ctx_set_decode_path": (_c_int, [_vp, _c_int]),
    "tq_quantize_kv": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _vp]),
    "tq_decode_workspace_bytes": (_c_size, [_vp, _c_int, _c_int, _c_int, _c_int]),
    "tq_attn_decode": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp, _vp,
                                _c_size, _vp]),
    "tq_attn_decode_noalloc": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp, _vp]),
    "tq_dequantize_kv": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp, _vp]),
    "tq_ip_topk_workspace_bytes": (_c_size, [_vp, _c_int, _c_int, _c_int, _c_int]),
    "tq_ip_topk": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _c_size,
                            _vp]),
    "tq_ctx_set_sparse_v": (_c_int, [_vp, ctypes.c_float]),
    "tq_paged_pool_bytes": (_c_size, [_vp, _c_int, _c_int]),
    "tq_quantize_kv_paged": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _c_int, _vp, _c_int, _vp]),
    "tq_attn_decode_paged": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _c_int, _vp, _vp, _vp,
                                      _vp, _c_size, _vp]),
    "tq_dequantize_kv_paged": (_c_int, [_vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp,
                                        _vp]),
    "tq_ip_topk_paged": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _c_int, _vp, _c_int, _vp,
                                  _vp, _vp, _c_size, _vp]),
    "tq_quantize_kv_strided": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(ctypes.c_int64), _c_int, _c_int, _c_int, _vp,
                                        _vp, _c_int, _vp]),
    "tq_quantize_kv_paged_strided": (_c_int, [_vp, _vp, _vp, ctypes.POINTER(ctypes.c_int64), _c_int, _c_int, _c_int,
                                              _vp, _vp, _c_int, _vp, _c_int, _vp]),
    "tq_selftest_bounded_wait": (_c_int, [_vp, _vp]),
    "tq_get_device_status": (_c_int, [_vp, _vp]),
    "tq_status_string": (ctypes.c_char_p, [_c_int]),
}


class TQError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")


def header_functions():
    """Names of the functions ``include/tq.h`` declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_\w+)\s*\(", text)))


def lib():
    """Loads libtq.so once (building it in-tree with nvcc first if it is missing or older
    than its sources).  Raises if that fails."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            if not _build.up_to_date():
                _build.build()
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status):
    return lib().tq_status_string(int(status)).decode()


def _check(fn, rc):
    if rc != TQ_OK:
        raise TQError(fn, rc)


def _ptr(t):
    """Device (or host) address of a tensor, or None."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---- host-only set-up ------------------------------------------------------------------

def tq_make_codebook(d, levels):
    """(centroids [levels], boundaries [levels-1]) as lists of floats (fp64)."""
    c = (ctypes.c_double * levels)()
    t = (ctypes.c_double * max(levels - 1, 1))()
    _check("tq_make_codebook", lib().tq_make_codebook(d, levels, c, t))
    return list(c), list(t)[:levels - 1]


def tq_make_rotation(d, seed):
    """Pi as a flat row-major list of d*d floats."""
    buf = (ctypes.c_double * (d * d))()
    _check("tq_make_rotation", lib().tq_make_rotation(d, ctypes.c_uint64(seed), buf))
    return list(buf)


def tq_make_projection(m, d, seed):
    """S as a flat row-major list of m*d floats."""
    buf = (ctypes.c_double * (m * d))()
    _check("tq_make_projection", lib().tq_make_projection(m, d, ctypes.c_uint64(seed), buf))
    return list(buf)


# ---- raw C-ABI wrappers (pointers are ints or ctypes values) -------------------------------

def tq_ctx_create(d, bits, m, seed, device):
    out = ctypes.c_void_p()
    _check("tq_ctx_create", lib().tq_ctx_create(d, bits, m, ctypes.c_uint64(seed), device, ctypes.byref(out)))
    return out


def tq_ctx_create_kv(d, key_bits, value_bits, qjl, seed, device):
    out = ctypes.c_void_p()
    _check("tq_ctx_create_kv", lib().tq_ctx_create_kv(d, key_bits, value_bits, 1 if qjl else 0, ctypes.c_uint64(seed),
                                                      device, ctypes.byref(out)))
    return out


def tq_ctx_destroy(ctx):
    lib().tq_ctx_destroy(ctx)


def tq_page_bytes(ctx):
    return lib().tq_page_bytes(ctx)


def tq_cache_bytes(ctx, batch, kv_heads, max_tokens):
    return lib().tq_cache_bytes(ctx, batch, kv_heads, max_tokens)


def tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens):
    return lib().tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens)


def tq_quantize_kv(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, stream):
    return lib().tq_quantize_kv(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, stream)


def tq_attn_decode(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                   workspace, workspace_bytes, stream):
    return lib().tq_attn_decode(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out,
                                logits_out, workspace, workspace_bytes, stream)


def tq_attn_decode_noalloc(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out, stream):
    return lib().tq_attn_decode_noalloc(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out,
                                        logits_out, stream)


def tq_get_device_status(ctx, stream):
    return lib().tq_get_device_status(ctx, stream)


def tq_status_string(status):
    return status_string(status)


def tq_ctx_get_constants(ctx, d, bits, m):
    """dict(pi, s, ck, tk, cv, tv) of flat fp64 lists (the context's host copies)."""
    lk, lv = 2 ** (bits - 1), 2 ** bits
    bufs = dict(pi=(ctypes.c_double * (d * d))(), s=(ctypes.c_double * (m * d))(),
                ck=(ctypes.c_double * lk)(), tk=(ctypes.c_double * (lk - 1))(),
                cv=(ctypes.c_double * lv)(), tv=(ctypes.c_double * (lv - 1))())
    _check("tq_ctx_get_constants", lib().tq_ctx_get_constants(ctx, bufs["pi"], bufs["s"], bufs["ck"], bufs["tk"],
                                                              bufs["cv"], bufs["tv"]))
    return {k: list(v) for k, v in bufs.items()}


# ---- tensor-level convenience (still only marshalling) --------------------------------------

class Context:
    """One (d, bits, m, seed) context on one CUDA device; wraps the C-ABI calls for torch
    tensors.  Every method is asynchronous on the given (or current) stream.  With key_bits
    (and value_bits, qjl) the context has separate key and value widths (format version 2,
    tq_ctx_create_kv); bits is then ignored."""

    def __init__(self, d, bits=None, m=None, seed=0, device=0, decode_path="auto", key_bits=None,
                 value_bits=None, qjl=True):
        self.d, self.seed, self.device = d, seed, device
        if key_bits is not None:
            self.key_bits, self.value_bits, self.qjl = key_bits, value_bits, bool(qjl)
            self.bits, self.m = None, d if qjl else 0
            self._ctx = tq_ctx_create_kv(d, key_bits, value_bits, qjl, seed, device)
        else:
            self.bits, self.m = bits, d if m is None else m
            self._ctx = tq_ctx_create(d, bits, self.m, seed, device)
        if decode_path != "auto":
            self.set_decode_path(decode_path)

    def set_decode_path(self, path):
        """'auto', 'simt', 'mma', 'tc' or 'tc4' (TQ_DECODE_*); query workspace sizes afterwards."""
        code = DECODE_PATHS[path] if isinstance(path, str) else int(path)
        _check("tq_ctx_set_decode_path", lib().tq_ctx_set_decode_path(self._ctx, code))
        self.decode_path = path

    def set_sparse_v(self, threshold):
        """Sparse V: positions with p_t = exp(l_t - running max) below threshold add no value
        (0 = dense attention, the default)."""
        _check("tq_ctx_set_sparse_v", lib().tq_ctx_set_sparse_v(self._ctx, float(threshold)))
        self.sparse_v = float(threshold)

    def close(self):
        if self._ctx:
            tq_ctx_destroy(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._ctx

    @property
    def page_bytes(self):
        return tq_page_bytes(self._ctx)

    def cache_bytes(self, batch, kv_heads, max_tokens):
        return tq_cache_bytes(self._ctx, batch, kv_heads, max_tokens)

    def workspace_bytes(self, batch, q_heads, kv_heads, max_tokens):
        return tq_decode_workspace_bytes(self._ctx, batch, q_heads, kv_heads, max_tokens)

    def alloc_cache(self, batch, kv_heads, max_tokens):
        import torch
        n = self.cache_bytes(batch, kv_heads, max_tokens)
        if n == 0:
            raise TQError("tq_cache_bytes", TQ_EINVAL)
        return torch.empty(n, dtype=torch.uint8, device=f"cuda:{self.device}")

    def alloc_workspace(self, batch, q_heads, kv_heads, max_tokens):
        import torch
        n = self.workspace_bytes(batch, q_heads, kv_heads, max_tokens)
        if n == 0:
            raise TQError("tq_decode_workspace_bytes", TQ_EINVAL)
        return torch.empty(n, dtype=torch.uint8, device=f"cuda:{self.device}")

    def quantize_kv(self, k, v, start_pos, cache, max_tokens, stream=None):
        """k, v: bf16 [B, Hkv, n_tokens, d] contiguous; start_pos: int32 [B] on the device."""
        B, H, N, d = k.shape
        rc = tq_quantize_kv(self._ctx, _ptr(k), _ptr(v), B, H, N, _ptr(start_pos), _ptr(cache), max_tokens,
                            _stream_handle(stream))
        _check("tq_quantize_kv", rc)

    def dequantize_kv(self, cache, start_pos, batch, kv_heads, n_tokens, max_tokens, k_out=None, v_out=None,
                      stream=None):
        """Reconstructed keys / values (fp32 [B, Hkv, n_tokens, d]) of the slots from start_pos[b]."""
        rc = lib().tq_dequantize_kv(self._ctx, _ptr(cache), batch, kv_heads, max_tokens, _ptr(start_pos), n_tokens,
                                    _ptr(k_out), _ptr(v_out), _stream_handle(stream))
        _check("tq_dequantize_kv", rc)

    def attn_decode(self, q, cache, seq_lens, kv_heads, max_tokens, out, workspace, logits=None, stream=None):
        """q, out: fp32 [B, Hq, d]; seq_lens: int32 [B] on the device; logits: None or
        fp32 [B, Hq, max_tokens]."""
        B, Hq, d = q.shape
        rc = tq_attn_decode(self._ctx, _ptr(q), B, Hq, kv_heads, _ptr(cache), _ptr(seq_lens), max_tokens,
                            _ptr(out), _ptr(logits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream_handle(stream))
        _check("tq_attn_decode", rc)

    @staticmethod
    def _kv_strides(k, v):
        """int64[6] element strides (batch, kv head, token) of k and v, viewed as [B, H, T, d]
        with unit stride in d (a permuted view of a [B, T, H, d] projection output is fine)."""
        if k.shape != v.shape or k.stride(3) != 1 or v.stride(3) != 1:
            raise TQError("tq_quantize_kv_strided", TQ_EINVAL)
        st = (ctypes.c_int64 * 6)(*(k.stride()[:3] + v.stride()[:3]))
        return st

    def quantize_kv_strided(self, k, v, start_pos, cache, max_tokens, stream=None):
        """quantize_kv for k, v of logical shape [B, Hkv, n_tokens, d] with any strides (unit in d)."""
        B, H, N, d = k.shape
        rc = lib().tq_quantize_kv_strided(self._ctx, _ptr(k), _ptr(v), self._kv_strides(k, v), B, H, N,
                                          _ptr(start_pos), _ptr(cache), max_tokens, _stream_handle(stream))
        _check("tq_quantize_kv_strided", rc)

    def quantize_kv_paged_strided(self, k, v, start_pos, pool, n_blocks, block_table, stream=None):
        B, H, N, d = k.shape
        rc = lib().tq_quantize_kv_paged_strided(self._ctx, _ptr(k), _ptr(v), self._kv_strides(k, v), B, H, N,
                                                _ptr(start_pos), _ptr(pool), n_blocks, _ptr(block_table),
                                                block_table.shape[1], _stream_handle(stream))
        _check("tq_quantize_kv_paged_strided", rc)

    # ---- paged (block-table) cache: pool of blocks, each the kv_heads pages of 128 slots ----
    def alloc_pool(self, kv_heads, n_blocks):
        import torch
        n = lib().tq_paged_pool_bytes(self._ctx, kv_heads, n_blocks)
        if n == 0:
            raise TQError("tq_paged_pool_bytes", TQ_EINVAL)
        return torch.empty(n, dtype=torch.uint8, device=f"cuda:{self.device}")

    def quantize_kv_paged(self, k, v, start_pos, pool, n_blocks, block_table, stream=None):
        """k, v: bf16 [B, Hkv, n_tokens, d]; block_table: int32 [B, max_blocks] on the device."""
        B, H, N, d = k.shape
        rc = lib().tq_quantize_kv_paged(self._ctx, _ptr(k), _ptr(v), B, H, N, _ptr(start_pos), _ptr(pool), n_blocks,
                                        _ptr(block_table), block_table.shape[1], _stream_handle(stream))
        _check("tq_quantize_kv_paged", rc)

    def attn_decode_paged(self, q, pool, n_blocks, block_table, seq_lens, kv_heads, out, workspace, logits=None,
                          stream=None):
        """As attn_decode, on a block pool; the workspace is that of max_tokens = 128 * max_blocks."""
        B, Hq, d = q.shape
        rc = lib().tq_attn_decode_paged(self._ctx, _ptr(q), B, Hq, kv_heads, _ptr(pool), n_blocks, _ptr(block_table),
                                        block_table.shape[1], _ptr(seq_lens), _ptr(out), _ptr(logits), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream_handle(stream))
        _check("tq_attn_decode_paged", rc)

    def dequantize_kv_paged(self, pool, n_blocks, block_table, start_pos, batch, kv_heads, n_tokens, k_out=None,
                            v_out=None, stream=None):
        rc = lib().tq_dequantize_kv_paged(self._ctx, _ptr(pool), n_blocks, _ptr(block_table), block_table.shape[1],
                                          batch, kv_heads, _ptr(start_pos), n_tokens, _ptr(k_out), _ptr(v_out),
                                          _stream_handle(stream))
        _check("tq_dequantize_kv_paged", rc)

    def ip_topk_paged(self, q, pool, n_blocks, block_table, seq_lens, kv_heads, k, out_idx=None, out_score=None,
                      workspace=None, stream=None):
        """ip_topk on a block pool (block_table int32 [B, max_blocks] on the device)."""
        import torch
        B, Hq, d = q.shape
        T = 128 * block_table.shape[1]
        if out_idx is None:
            out_idx = torch.empty(B, Hq, k, dtype=torch.int32, device=q.device)
        if out_score is None:
            out_score = torch.empty(B, Hq, k, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = self.alloc_topk_workspace(B, Hq, kv_heads, T)
        rc = lib().tq_ip_topk_paged(self._ctx, _ptr(q), B, Hq, kv_heads, _ptr(pool), n_blocks, _ptr(block_table),
                                    block_table.shape[1], _ptr(seq_lens), k, _ptr(out_idx), _ptr(out_score),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream))
        _check("tq_ip_topk_paged", rc)
        return out_idx, out_score

    def alloc_topk_workspace(self, batch, q_heads, kv_heads, max_tokens, device="cuda"):
        """Device scratch of tq_ip_topk (tq_ip_topk_workspace_bytes bytes)."""
        import torch
        n = lib().tq_ip_topk_workspace_bytes(self._ctx, batch, q_heads, kv_heads, max_tokens)
        if n == 0:
            raise TQError("tq_ip_topk_workspace_bytes", TQ_EINVAL)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def ip_topk(self, q, cache, seq_lens, kv_heads, max_tokens, k, out_idx=None, out_score=None, workspace=None,
                stream=None):
        """Compressed inner-product scan (tq_ip_topk): per query head the k slots with the largest
        estimated <q, k^_t>.  q: fp32 [B, Hq, d]; seq_lens: int32 [B] on the device.  Returns
        (out_idx int32 [B, Hq, k], out_score fp32 [B, Hq, k])."""
        import torch
        B, Hq, d = q.shape
        if out_idx is None:
            out_idx = torch.empty(B, Hq, k, dtype=torch.int32, device=q.device)
        if out_score is None:
            out_score = torch.empty(B, Hq, k, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = self.alloc_topk_workspace(B, Hq, kv_heads, max_tokens)
        rc = lib().tq_ip_topk(self._ctx, _ptr(q), B, Hq, kv_heads, _ptr(cache), _ptr(seq_lens), max_tokens, k,
                              _ptr(out_idx), _ptr(out_score), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream))
        _check("tq_ip_topk", rc)
        return out_idx, out_score

    def device_status(self, stream=None):
        """Synchronises the stream; returns (and clears) the sticky device status code."""
        return tq_get_device_status(self._ctx, _stream_handle(stream))

    def constants(self):
        return tq_ctx_get_constants(self._ctx, self.d, self.bits, self.m)
