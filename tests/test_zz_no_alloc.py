"""The allocation-free split-KV call against the workspace call, through the C ABI.

mslk_attn_split_kv_static runs the same split-KV path as mslk_attn_split_kv but keeps its
workspace in a fixed array inside the library, for callers that cannot allocate device
memory when they call.  This file is collected after the other test files, so a run that
stops at the first failure has run everything else first; it also passes on its own.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

import attention_fmha_fwd_gb300 as fa
from attention_fmha_fwd_gb300 import _capi, build, inputs
from tests.gpu_util import compare


def test_static_workspace_limit_is_enforced_before_launch():
    """A problem whose workspace exceeds the fixed array is refused with a reason before
    anything is launched (no GPU needed)."""
    build.build()
    lib = _capi.load()
    a = _capi.AttnArgs()
    a.q = a.k = a.v = a.out = a.lse = 0x10000  # never dereferenced: the size check comes first
    a.B, a.M, a.Mkv, a.H, a.Hkv, a.K, a.Kv = 8, 1024, 8192, 16, 0, 128, 128
    a.sq = a.so = _capi.Strides(1024 * 16 * 128, 16 * 128, 128)
    a.sk = a.sv = _capi.Strides(8192 * 16 * 128, 16 * 128, 128)
    # 64 chunks of fp32 [8, 1024, 16, 128] outputs: 4 GiB, far beyond the fixed array
    st = lib.mslk_attn_split_kv_static(ctypes.byref(a), 64, None)
    assert st == _capi.MSLK_ERR_UNSUPPORTED
    why = lib.mslk_last_error().decode()
    assert "fixed" in why and str(_capi.SPLIT_KV_STATIC_BYTES) in why


@pytest.mark.gpu
def test_static_split_kv_matches_workspace_call_twice():
    """Two calls in a row (different problems, so the second finds the first's data in the
    array): each equals the workspace call within the parity tolerances, and neither
    allocates device memory."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    cases = [(1, 128, 1024, 16, 128, 8, "none", {}),           # the split-KV workload
             (2, 200, 1500, 4, 64, 5, "causal_bottom_right", {})]
    for B, M, Mkv, H, D, n, mask, kw in cases:
        q, k, v = (t.cuda() for t in inputs.qkv(B, M, Mkv, H, D, seed=60 + n))
        ref_out, ref_lse = fa.attn_split_kv(q, k, v, n_chunks=n, mask=mask, **kw)
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        torch.cuda.synchronize()
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        fa.attn_split_kv_static(q, k, v, n_chunks=n, mask=mask, out=out, lse=lse, **kw)
        torch.cuda.synchronize()
        assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == before
        compare(out.double().cpu().numpy(), lse.double().cpu().numpy(),
                ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                f"static split B{B} M{M} Mkv{Mkv} n{n} {mask}")
    assert fa.device_status() == 0
