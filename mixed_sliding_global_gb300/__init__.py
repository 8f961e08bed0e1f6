"""Mixed sliding/global GQA attention over a device-resident KV cache, for NVIDIA GB300.

Python binding of the C ABI in ``include/gemma_attn.h`` (``libgemma_attn.so``). The functions
below carry the C names and only marshal arguments: sizes are read from tensor shapes,
pointers from ``data_ptr()``, and the stream from torch's current stream. Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
loading fails loudly when the library has not been built.
"""
from .binding import (  # noqa: F401
    GEMMA_SLIDING, GEMMA_GLOBAL, GEMMA_SLIDING_RING, GEMMA_BF16, GEMMA_FP32, GEMMA_OK,
    GEMMA_DEVERR_SEQ_LEN, GEMMA_DEVERR_WRITE_POS, GEMMA_DEVERR_TIMEOUT, GEMMA_DEVERR_N_REAL,
    GEMMA_DEVERR_PAGE,
    GemmaError, library, library_path, exported_symbols,
    gemma_kv_append, gemma_attn_decode, gemma_attn_decode_static, gemma_attn_prefill, gemma_attn_softcap,
    gemma_kv_append_bucket, gemma_attn_prefill_bucket, gemma_attn_decode_append,
    gemma_kv_append_ring, gemma_kv_append_paged, gemma_attn_paged, gemma_attn_workspace_size_paged,
    gemma_attn_workspace_size, gemma_logit_softcap_argmax, gemma_logit_workspace_size,
    gemma_status_string, gemma_abi_version,
)
