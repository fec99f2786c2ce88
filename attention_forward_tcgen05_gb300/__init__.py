"""GB300 (sm_103a) attention-forward engine: exact SDPA with online softmax.

Prefill FMHA on tcgen05 tensor cores (TMA-fed, TMEM accumulators) and a GQA
split-KV decode with an LSE-weighted merge, behind the C ABI of
``include/attn.h``.  ``libattn.so`` is built in-tree by ``build.build()``.
"""
from ._binding import (  # noqa: F401
    ATTN_BF16, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_INPUT, ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_INVALID_ARG,
    ATTN_ERR_SCRATCH_TOO_SMALL, ATTN_ERR_UNSUPPORTED, ATTN_F32, ATTN_OK, LIB_PATH, AttnError,
    attn_debug_wait_timeout, attn_decode, attn_decode_noalloc, attn_decode_noalloc_scratch_bytes,
    attn_decode_packed, attn_decode_split, attn_decode_split_packed, attn_merge, attn_prefill_fwd,
    attn_prefill_packed, attn_prefill_schedule, attn_prefill_varlen, attn_prefill_varlen_window,
    attn_prefill_window, attn_strerror, attn_sync_check, attn_version, decode, decode_counters,
    decode_packed, decode_split, decode_split_packed, load, merge, prefill, prefill_schedule,
    prefill_varlen, prefill_window, sync_check)
