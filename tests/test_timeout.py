"""Bounded waits: a wait nobody signals ends with an error status, not a hang."""
import ctypes

import pytest
import torch

import attention_forward_tcgen05_gb300 as attn

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_context_survives():
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert attn.attn_sync_check(s) == attn.ATTN_OK
    assert attn.attn_debug_wait_timeout(2_000_000, s) == attn.ATTN_OK  # 2 ms limit
    assert attn.attn_sync_check(s) == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_sync_check(s) == attn.ATTN_OK  # the error word was cleared
    # the context is still usable
    q = torch.randn(1, 130, 2, 64, device="cuda").to(torch.bfloat16)
    o, lse = attn.prefill(q, q, q, causal=True)
    assert attn.attn_sync_check(s) == attn.ATTN_OK
    assert torch.isfinite(o.float()).all()
