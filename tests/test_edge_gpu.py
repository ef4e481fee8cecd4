"""Numerical and shape edge cases on both kernels, vs the fp64 oracle through the C ABI.

* large logits (scale x 30: scores hundreds apart), so the lazy rescale and the empty
  -inf handling work at the extremes of fp32 exponents;
* a key late in the row that dominates it (the running max jumps after many tiles);
* many key tiles per row (accumulation over 512 tiles, sampled rows);
* unit counts that do not divide the SM count, and many heads on the decode path.
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

KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL}


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


def _run(q, k, v, scale, mask, policy=0):
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=scale)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("M,Mkv,mask,policy", [
    (300, 900, "none", 0), (300, 300, "causal", 0), (4, 3000, "none", 0), (4, 3000, "none", 1)])
def test_large_logits(M, Mkv, mask, policy):
    """scale 30/sqrt(D): logits span hundreds; softmax is near one-hot per row."""
    q, k, v = inputs.qkv(1, M, Mkv, 2, 128, seed=M + Mkv)
    s = 30.0 / 128 ** 0.5
    out, lse = _run(q, k, v, s, mask, policy)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask])
    compare(out, lse, ro, rl, f"large logits M{M} Mkv{Mkv} {mask} policy{policy}")


@pytest.mark.parametrize("M,policy", [(256, 0), (2, 0), (2, 1)])
def test_late_dominant_key(M, policy):
    """Key Mkv - 5 has a large dot product with every query: the running max jumps by far
    more than the lazy threshold in the last tile, after many tiles of small scores."""
    Mkv, H, D = 4000, 2, 128
    q, k, v = inputs.qkv(1, M, Mkv, H, D, seed=41)
    k = k.clone()
    qm = q.float().mean(dim=1, keepdim=True)            # [1, 1, H, D]
    k[:, Mkv - 5] = (qm[:, 0] * 40.0).to(torch.bfloat16)  # aligned with the average query
    s = D ** -0.5
    out, lse = _run(q, k, v, s, "none", policy)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out, lse, ro, rl, f"late dominant key M{M} policy{policy}")


def test_many_key_tiles_sampled():
    """256 queries against 65536 keys (512 key tiles per row), rows sampled for the oracle."""
    M, Mkv, H, D = 256, 65536, 2, 128
    q, k, v = inputs.qkv(1, M, Mkv, H, D, seed=8)
    s = D ** -0.5
    out, lse = _run(q, k, v, s, "causal")  # top-left causal: row i sees keys 0..i
    out2, lse2 = fa.attn_fwd(*to_dev(q, k, v), mask="none", scale=s)
    out2, lse2 = out2.double().cpu().numpy(), lse2.double().cpu().numpy()
    rows = [0, 1, 77, 128, 255]
    qs = q[:, rows]
    ro, rl = oracle.attention(f32(qs), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out2[:, rows], lse2[:, :, rows], ro, rl, "65536 keys, sampled rows")
    # causal: row i against its own prefix
    for i in (0, 77, 255):
        ro, rl = oracle.attention(f32(q[:, i:i + 1]), f32(k[:, :i + 1]), f32(v[:, :i + 1]), s,
                                  oracle.MASK_NONE)
        compare(out[:, i:i + 1], lse[:, :, i:i + 1], ro, rl, f"causal row {i}")


@pytest.mark.parametrize("B,M,Mkv,H,D,mask", [
    (3, 300, 300, 40, 64, "causal"),     # 3 x 40 x 2 = 240 units on 152 SMs
    (5, 1, 1000, 96, 128, "none"),       # 480 decode CTAs
    (1, 7, 513, 128, 64, "causal"),      # 128 heads, 7 rows
])
def test_odd_unit_counts(B, M, Mkv, H, D, mask):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=B * H + M)
    s = D ** -0.5
    out, lse = _run(q, k, v, s, mask)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask])
    compare(out, lse, ro, rl, f"B{B} M{M} Mkv{Mkv} H{H} D{D} {mask}")


@pytest.mark.parametrize("M,policy", [(4, 0), (4, 2), (8, 0), (2, 0)])
def test_few_rows_many_heads_dispatch(M, policy):
    """Few query rows over 16 x 8 (batch, head) units: the automatic choice sends 2+ rows to
    the tensor cores (policy 0), policy 2 keeps the CUDA-core kernel; both match the oracle."""
    B, Mkv, H, D = 16, 3000, 8, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=M + 100)
    s = D ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="causal", scale=s, bottom_right=True)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_CAUSAL, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"M{M} policy{policy}")
