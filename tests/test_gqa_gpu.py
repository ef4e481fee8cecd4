"""Grouped-query attention (Hkv K/V heads for H query heads): CUDA path vs the fp64 oracle.

Query head h reads K/V head h // (H / Hkv) (the pages' BMGHK layout flattened group-major).
Few query rows fold a group's query heads into one block of rows (each K/V head streamed
once); the tensor-core path maps heads per unit.  All calls go through the C ABI
(mslk_attn with Hkv set).
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

KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL,
        "blockdiag": oracle.MASK_BLOCKDIAG, "blockdiag_causal": oracle.MASK_BLOCKDIAG_CAUSAL}


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


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def _np(t):
    return t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


@pytest.mark.parametrize("B,M,Mkv,H,Hkv,D,mask,br,wl,policy", [
    (2, 1, 3000, 8, 2, 128, "causal", True, None, 0),     # decode, 4 heads folded per K/V head
    (1, 2, 2500, 8, 2, 128, "causal", True, None, 0),     # 2 positions x 4 heads = 8 rows
    (1, 3, 2000, 8, 2, 64, "causal", True, 100, 0),       # 3 positions: 2 heads folded
    (2, 4, 1500, 6, 3, 128, "none", False, None, 0),      # group 2, 4 positions: 2 heads folded
    (1, 1, 5000, 16, 1, 128, "none", False, None, 0),     # one K/V head for 16 query heads (fold 8)
    (1, 300, 700, 8, 2, 128, "causal", True, None, 0),    # tensor cores
    (2, 260, 260, 6, 2, 64, "causal", False, 50, 0),
    (1, 4, 900, 8, 4, 128, "causal", True, None, 1),      # few rows forced onto the tensor cores
])
def test_gqa_dense(B, M, Mkv, H, Hkv, D, mask, br, wl, policy):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, Hkv=Hkv, seed=M + H + Hkv)
    s = D ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=br, window_left=wl)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=br, window_left=wl)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"gqa B{B} M{M} Mkv{Mkv} H{H}/{Hkv} D{D} {mask} policy{policy}")


@pytest.mark.parametrize("lq", [[1, 1, 1], [2, 1, 2], [100, 7, 300]])
def test_gqa_varlen(lq):
    lk = [900, 64, 1300]
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q, k, v = inputs.qkv(1, sum(lq), sum(lk), 8, 128, Hkv=2, seed=sum(lq))
    s = 128 ** -0.5
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", scale=s, cu_seqlens_q=_i32(cu_q),
                           cu_seqlens_k=_i32(cu_k), max_seqlen_q=max(lq), max_seqlen_k=max(lk),
                           bottom_right=True)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k,
                              bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"gqa varlen {lq}")


def test_gqa_paged_decode():
    lq, lk, ps, H, Hkv = [1, 1, 2], [700, 3001, 129], 64, 8, 2
    table, n_pages, _ = inputs.page_table(lk, ps, spare_pages=2, seed=4)
    q, k, v = inputs.qkv(1, sum(lq), n_pages * ps, H, 128, Hkv=Hkv, seed=4)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd_lanes(q.cuda(), k.cuda().view(n_pages, ps, Hkv, 128),
                                 v.cuda().view(n_pages, ps, Hkv, 128), seqlen_k=_i32(lk),
                                 cu_seqlens_q=_i32(inputs.cu_seqlens(lq)), max_seqlen_q=max(lq),
                                 max_seqlen_k=max(lk), block_table=table.cuda(), page_size=ps,
                                 bottom_right=True)
    ro, rl = oracle.attention_lanes(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL,
                                    inputs.cu_seqlens(lq), lk, block_table=table.numpy(),
                                    page_size=ps, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "gqa paged decode")


@pytest.mark.parametrize("M", [1, 200])
def test_gqa_split_kv(M):
    q, k, v = inputs.qkv(2, M, 2048, 8, 128, Hkv=2, seed=M)
    s = 128 ** -0.5
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in inputs.equal_chunks(2048, 4):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=s, kv_offset=a)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"gqa split-KV M{M}")


def test_gqa_fp8_decode():
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(2, 1, 4000, 8, 128, Hkv=2, seed=3)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(),
                               mask="causal", scale=s, bottom_right=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), s,
                                  oracle.MASK_CAUSAL, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "gqa fp8 decode")


def test_gqa_equals_expanded_on_tensor_cores():
    """Grouped heads give the same bits as the same K/V repeated per query head (the tensor
    cores process each query head's unit the same way in both)."""
    q, k, v = inputs.qkv(1, 400, 400, 8, 128, Hkv=2, seed=17)
    qd, kd, vd = to_dev(q, k, v)
    a = fa.attn_fwd(qd, kd, vd, mask="causal")
    b = fa.attn_fwd(qd, kd.repeat_interleave(4, dim=2), vd.repeat_interleave(4, dim=2), mask="causal")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ folded heads on the tensor cores
# One query position per batch / sequence, group > 1, and >= 64 (batch, K/V head) units
# (or the tensor-core policy): the group's query heads become the rows of one unit.

@pytest.mark.parametrize("B,Mkv,H,Hkv,D,mask,br,wl,policy", [
    (16, 3000, 32, 4, 128, "causal", True, None, 0),     # 64 units, bottom-right causal
    (8, 2500, 64, 8, 64, "causal", True, 200, 0),        # window relative to the last key
    (16, 700, 16, 4, 128, "causal", False, None, 0),     # top-left: the query sees key 0 only
    (2, 2000, 24, 2, 128, "none", False, None, 1),       # few units, forced onto the tensor cores
    (64, 300, 16, 1, 128, "none", False, None, 0),       # one K/V head for 16 query heads
])
def test_folded_heads_dense(B, Mkv, H, Hkv, D, mask, br, wl, policy):
    q, k, v = inputs.qkv(B, 1, Mkv, H, D, Hkv=Hkv, seed=B + Mkv + H)
    s = D ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=br, window_left=wl)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=br, window_left=wl)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"folded B{B} Mkv{Mkv} H{H}/{Hkv} D{D} {mask} br{br} wl{wl}")


def test_folded_heads_varlen_and_paged():
    """70 packed sequences with one query each (some with none), 2 K/V heads of 4 query heads."""
    n = 70
    g = torch.Generator().manual_seed(12)
    lq = [0 if i % 9 == 4 else 1 for i in range(n)]
    lk = torch.randint(1, 1500, (n,), generator=g).tolist()
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q, k, v = inputs.qkv(1, sum(lq), sum(lk), 8, 128, Hkv=2, seed=12)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", scale=s, cu_seqlens_q=_i32(cu_q),
                           cu_seqlens_k=_i32(cu_k), max_seqlen_q=1, max_seqlen_k=max(lk),
                           bottom_right=True)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k,
                              bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "folded varlen")
    # the same lanes paged (128-key pages)
    ps = 128
    table, n_pages, _ = inputs.page_table(lk, ps, spare_pages=1, seed=12)
    rows = np.concatenate([oracle.lane_rows(i, lk, block_table=table.numpy(), page_size=ps) for i in range(n)])
    kp = torch.zeros((1, n_pages * ps, 2, 128), dtype=torch.bfloat16)
    vp = torch.zeros((1, n_pages * ps, 2, 128), dtype=torch.bfloat16)
    kp[0, torch.from_numpy(rows)] = k[0]
    vp[0, torch.from_numpy(rows)] = v[0]
    out, lse = fa.attn_fwd_lanes(q.cuda(), kp.cuda().view(n_pages, ps, 2, 128),
                                 vp.cuda().view(n_pages, ps, 2, 128), seqlen_k=_i32(lk),
                                 cu_seqlens_q=_i32(cu_q), max_seqlen_q=1, max_seqlen_k=max(lk),
                                 block_table=table.cuda(), page_size=ps, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "folded paged")


def test_folded_heads_partial_merge():
    q, k, v = inputs.qkv(32, 1, 2048, 16, 128, Hkv=2, seed=21)
    s = 128 ** -0.5
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in inputs.equal_chunks(2048, 3):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=s, mask="causal", kv_offset=a - 2047)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_CAUSAL, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "folded split-KV")


def test_folded_heads_fp8():
    """E4M3 with per-head descales: every folded row has its own query descale."""
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(16, 1, 2500, 16, 128, Hkv=4, seed=5)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(),
                               mask="causal", scale=s, bottom_right=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), s,
                                  oracle.MASK_CAUSAL, bottom_right=True)
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.abs(lse - rl).max() <= 1e-3
    # E4M3 probabilities on the tensor cores: |d out| <= 2^-4 sum p|v| / sum p (+ output rounding)
    from tests.test_fp8_gpu import _deq, _p_rounding_check
    _p_rounding_check(out, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), s, "causal",
                      "folded fp8", br=True)
