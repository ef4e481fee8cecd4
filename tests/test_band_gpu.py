"""Bottom-right alignment and local windows: CUDA path vs the fp64 oracle, through the C ABI.

Masks of "Attention - Biases & masks" (LowerTriangularFromBottomRightMask, the local
attention masks, the block-diagonal bottom-right and local variants), in the reading the
oracle documents: query i pairs with key i + (bottom_right ? Lk - Lq : 0); windows keep
window_left keys before and window_right keys after the paired key.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fmha_fwd_gb300 as fa
import oracle
from attention_fmha_fwd_gb300 import inputs
from tests.gpu_util import compare, f32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_fmha_fwd_gb300 import build
    build.build()
    fa.set_path_policy(0)
    yield
    fa.set_path_policy(0)
    assert fa.device_status() == 0


KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL}


def _dense(B, M, Mkv, H, D, mask, br=False, wl=None, wr=None, seed=0, policy=0):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=seed)
    s = 1 / D ** 0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=br,
                               window_left=wl, window_right=wr)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=br,
                              window_left=wl, window_right=wr)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"B{B} M{M} Mkv{Mkv} H{H} D{D} {mask} br{br} wl{wl} wr{wr} policy{policy}")


@pytest.mark.parametrize("B,M,Mkv,H,D,mask,br,wl,wr", [
    (1, 300, 700, 2, 128, "causal", True, None, None),     # bottom-right causal, Mkv > M
    (2, 500, 200, 2, 64, "causal", True, None, None),      # M > Mkv: leading rows see nothing
    (1, 777, 777, 2, 128, "causal", False, 100, None),     # causal window, tiles skipped
    (1, 256, 1000, 2, 128, "causal", True, 63, None),      # bottom-right causal window
    (1, 600, 650, 2, 64, "none", True, 130, 70),           # two-sided local window
    (1, 300, 300, 2, 128, "none", False, 0, 0),            # one key per row
    (1, 400, 900, 3, 128, "none", False, None, 40),        # right edge only
    (1, 1100, 1100, 2, 128, "causal", False, 300, None),   # several units, window < unit
])
def test_band_tensor_core(B, M, Mkv, H, D, mask, br, wl, wr):
    _dense(B, M, Mkv, H, D, mask, br, wl, wr, seed=M + Mkv)


@pytest.mark.parametrize("M,Mkv,mask,br,wl,wr", [
    (1, 3000, "causal", True, None, None),
    (5, 3000, "causal", True, 200, None),
    (8, 2500, "none", True, 100, 3),
    (3, 5000, "causal", False, None, None),    # top-left: only keys 0..2
    (7, 40000, "causal", True, 20000, None),   # long window: cluster split of the band
])
def test_band_decode_and_both_paths(M, Mkv, mask, br, wl, wr):
    _dense(2, M, Mkv, 2, 128, mask, br, wl, wr, seed=M, policy=2)   # CUDA-core kernel
    _dense(2, M, Mkv, 2, 128, mask, br, wl, wr, seed=M, policy=1)   # tensor-core kernel


@pytest.mark.parametrize("br,wl", [(True, None), (False, 64), (True, 100)])
def test_band_blockdiag(br, wl):
    """Packed sequences with unequal query and key lengths per sequence."""
    lq, lk = [100, 300, 50, 260], [200, 300, 400, 129]
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q, k, v = inputs.qkv(1, sum(lq), sum(lk), 2, 128, seed=9)
    s = 1 / 128 ** 0.5
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", scale=s, cu_seqlens_q=cq,
                           cu_seqlens_k=ck, max_seqlen_q=max(lq), max_seqlen_k=max(lk),
                           bottom_right=br, window_left=wl)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k,
                              bottom_right=br, window_left=wl)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"blockdiag br{br} wl{wl}")


def test_bottom_right_mask_kinds():
    """The shorthand kinds 4/5 equal causal + bottom_right."""
    q, k, v = inputs.qkv(1, 200, 450, 2, 64, seed=4)
    a = fa.attn_fwd(*to_dev(q, k, v), mask="causal_bottom_right")
    b = fa.attn_fwd(*to_dev(q, k, v), mask="causal", bottom_right=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    lq, lk = [70, 130], [150, 200]
    cq = torch.tensor(inputs.cu_seqlens(lq), dtype=torch.int32, device="cuda")
    ck = torch.tensor(inputs.cu_seqlens(lk), dtype=torch.int32, device="cuda")
    q, k, v = inputs.qkv(1, 200, 350, 2, 64, seed=5)
    kw = dict(cu_seqlens_q=cq, cu_seqlens_k=ck, max_seqlen_q=130, max_seqlen_k=200)
    a = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal_bottom_right", **kw)
    b = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", bottom_right=True, **kw)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("M", [4, 640])
def test_windowed_split_kv(M):
    """A causal window over chunks: windowed partials (kv_offset per chunk) merged equal the
    windowed forward of the oracle."""
    q, k, v = inputs.qkv(1, M, 1024, 2, 128, seed=12)
    s = 1 / 128 ** 0.5
    off = 1024 - M  # bottom-right alignment folded into kv_offset
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in ((0, 300), (300, 700), (700, 1024)):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], mask="causal", scale=s,
                                kv_offset=a - off, window_left=256)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_CAUSAL, bottom_right=True,
                              window_left=256)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"windowed split M{M}")
