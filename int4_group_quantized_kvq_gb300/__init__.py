"""INT4 group-quantized paged KV cache for NVIDIA GB300 (sm_103a).

The compute lives in ``libkvq.so`` (hand-written CUDA kernels behind the C ABI of
``include/kvq.h``); this package is its ctypes binding.  PyTorch is used only for
device memory and streams.

    from int4_group_quantized_kvq_gb300 import config, kvq_pool_bytes, kvq_quantize_append, ...
"""
from .binding import (  # noqa: F401
    ABI_SYMBOLS,
    KVQ_EINVAL,
    KVQ_ECUDA,
    KVQ_EUNSUPPORTED,
    KVQ_EWORKSPACE,
    KVQ_FLAG_BAD_PAGE,
    KVQ_FLAG_BAD_POSITION,
    KVQ_FLAG_WAIT_TIMEOUT,
    KVQ_OK,
    CacheConfig,
    KvqError,
    config,
    kvq_block_bytes,
    kvq_decode_attention,
    kvq_decode_attention_noalloc,
    kvq_decode_attention_window,
    kvq_decode_step,
    kvq_decode_step_window,
    kvq_decode_workspace_bytes,
    kvq_dequantize_to_fp16_pool,
    kvq_fp16_append,
    kvq_fp16_decode_attention,
    kvq_fp16_decode_workspace_bytes,
    kvq_fp16_pool_bytes,
    kvq_int8_decode_attention,
    kvq_int8_decode_workspace_bytes,
    kvq_int8_pool_bytes,
    kvq_int8_quantize_append,
    kvq_mixed_decode_attention,
    kvq_mixed_decode_workspace_bytes,
    new_fp16_workspace,
    kvq_dequantize,
    kvq_last_error,
    kvq_pool_bytes,
    kvq_quantize_append,
    kvq_read_status,
    kvq_version,
    lib,
    new_workspace,
)
