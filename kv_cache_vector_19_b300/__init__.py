"""TurboQuant compressed KV cache for one B300 (sm_103a): online quantizer + decode attention.

The compute path is ``libtq.so`` (CUDA kernels behind the C ABI in ``include/tq.h``);
``binding`` is its ctypes shim and ``workloads`` draws seeded synthetic inputs.
"""
from .binding import (DECODE_PATHS, PAGE_TOKENS, TQ_DECODE_AUTO, TQ_DECODE_MMA, TQ_DECODE_SIMT, TQ_DECODE_TC,
                      TQ_EBOUNDS, TQ_ECUDA, TQ_EINVAL, TQ_ENOMEM, TQ_ENOTCONV, TQ_ESCRATCH, TQ_ETIMEOUT,
                      TQ_EUNSUPPORTED, TQ_OK, Context, TQError, lib, tq_attn_decode,
                      tq_attn_decode_noalloc, tq_cache_bytes, tq_ctx_create, tq_ctx_destroy, tq_ctx_get_constants,
                      tq_decode_workspace_bytes, tq_get_device_status, tq_make_codebook, tq_make_projection,
                      tq_make_rotation, tq_page_bytes, tq_quantize_kv, tq_status_string)
