"""Failure detection without a GPU fault: a bounded in-kernel wait that runs out ends the
kernel cleanly, the host reads MSLK_ERR_DEVICE_TIMEOUT, and the context stays usable."""

import pytest
import torch

import attention_fmha_fwd_gb300 as fa
from attention_fmha_fwd_gb300 import _capi, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert fa.device_status() == _capi.MSLK_OK
    fa.set_wait_timeout_ns(200_000_000)  # 0.2 s
    try:
        fa.diag_bounded_wait()          # waits on a barrier nothing completes
        assert fa.device_status() == _capi.MSLK_ERR_DEVICE_TIMEOUT
        assert "bounded wait" in fa.last_error()
        assert fa.device_status() == _capi.MSLK_OK  # the word was cleared
    finally:
        fa.set_wait_timeout_ns(2_000_000_000)
    # the device still computes
    q, k, v = inputs.qkv(1, 64, 64, 1, 64, seed=0)
    out, lse = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert fa.device_status() == _capi.MSLK_OK
