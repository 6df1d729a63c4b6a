"""Failure paths on the GPU without faulting it: a bounded wait that runs
out, and host validation that refuses bad arguments before any launch."""

import pytest
import torch

from exact_tiled_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_timeout_reported_and_context_survives(fa):
    assert fa.fa_device_status() == fa.FA_OK
    assert fa.fa_selftest_wait_timeout(50_000_000) == fa.FA_OK  # 50 ms
    assert fa.fa_device_status(clear=True) == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status() == fa.FA_OK
    q, k, v = W.dense_inputs(1, 130, 2, 64, 5, "cuda")
    o, lse = fa.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_invalid_arguments_rejected(fa):
    q, k, v = W.dense_inputs(1, 64, 2, 64, 6, "cuda")
    o = torch.empty_like(q)
    assert fa.fa_fwd(q, k, v, o, None, 1, 2, 2, 64, 80, 0.1, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd(q, k, v, o, None, 1, 2, 2, 64, 64, -1.0, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(q, k, v, o, None, 1, 2, 3, 64, 64, 0.1, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(q.data_ptr() + 2, k, v, o, None, 1, 2, 2, 64, 64, 0.1, 0) == fa.FA_ERR_INVALID
    assert fa.fa_device_status() == fa.FA_OK
